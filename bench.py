"""Benchmark of the Fathom decode step on GB300.

One step = one decode step over all layers of the workload: per layer, the
per-query-group plan, the gather of the planned plane runs (host-resident
regime), the scan + top-k and the exact sparse attention over the winners,
for every (sequence, KV head) unit of the layer.  The reported value is
microseconds per layer-step (whole job: time / (steps * layers * sessions));
the JSON line also carries the scanned-bytes rate, the roofline of the
dominant kernel, the end-to-end figure through the C ABI with host buffers,
the clocks seen and the CPU oracle baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload host_1m]
                    [--budget 48] [--impl fathom|reference] [--fixed]

Multi-GPU: one process per GPU (torchrun); every rank serves its own session
(its own seeded store), no data-path collective ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_plane_kv_gb300 import synth  # noqa: E402

METRIC = "decode-step µs/layer and scan GB/s (% of PCIe/HBM roofline) at 1M tokens"
CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if torch.cuda.is_available() and local < torch.cuda.device_count():
        torch.cuda.set_device(local)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The largest of the ranks' values (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(w: synth.Workload, rank: int) -> synth.Workload:
    """Every rank serves its own session: the same shapes with a rank-specific seed
    (rank 0 keeps the workload's own seed).  Units are never split across ranks."""
    return synth.shrink(w, seed=w.seed + 1000003 * rank) if rank else w


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling every 10 ms with timestamps; stop() keeps the samples that fall
    inside the timed region (host wall-clock window), or, when the region is shorter than
    the sampling period, the samples nearest to it."""

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self, wait_s=3.0):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "10"], stdout=self.fh, stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < wait_s and os.path.getsize(self.path) == 0:
                time.sleep(0.02)
        except Exception:
            self.proc = None

    @staticmethod
    def _epoch(ts):
        import datetime
        try:
            return datetime.datetime.strptime(ts.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self, device_index=0, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.03)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10 or not f[1].isdigit() or int(f[1]) != device_index:
                continue
            rows.append((self._epoch(f[0]), f[1:]))
        os.unlink(self.path)
        inside = rows
        how = "all samples"
        if window and rows and all(t is not None for t, _ in rows):
            a, b = window
            inside = [r for r in rows if a <= r[0] <= b]
            how = "inside the timed region"
            if not inside:   # region shorter than the sampling period: the nearest samples
                rows.sort(key=lambda r: min(abs(r[0] - a), abs(r[0] - b)))
                inside = rows[:2]
                how = "nearest to the timed region (shorter than the 10 ms period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for _, r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for _, r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, r in inside for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": how}


# ---------------------------------------------------------------- workload
class Setup:
    """Builds the store and rows of one session on this rank (untimed)."""

    def __init__(self, w: synth.Workload, budget: int, rank: int, steps_total: int, fixed: bool,
                 path: str = "fused", groups: int = 4, want_theta: bool = False):
        from bit_plane_kv_gb300 import binding as B
        self.B = B
        self.w, self.budget, self.fixed = w, budget, fixed
        # the decode step needs the depths and the run list; theta (the water level)
        # is a diagnostic, requested only with --plan-theta
        self.want_theta = want_theta
        w = rank_workload(w, rank)
        self.L, self.H = w.layers, w.units_per_layer()
        self.n, self.G, self.D, self.k = w.n, w.G, w.D, w.k
        self.nb = B.nblocks(self.n)
        self.host = w.regime == "host"
        self.shape = B.make_shape(self.H, self.n, self.D, self.G, self.k, w.n_sink, w.n_recent)
        dev = "cuda"
        L, H, n, D, nb = self.L, self.H, self.n, self.D, self.nb
        t0 = time.time()
        alloc = (lambda *s, dtype: torch.empty(*s, dtype=dtype, pin_memory=True)) if self.host else \
                (lambda *s, dtype: torch.empty(*s, dtype=dtype, device=dev))
        self.planes = alloc(L, H, D, 4, nb, dtype=torch.int64)
        self.scales = alloc(L, H, D, nb, dtype=torch.int16)
        self.krows = alloc(L, H, n, D, dtype=torch.bfloat16)
        self.vrows = alloc(L, H, n, D, dtype=torch.bfloat16)
        self.var = torch.empty(L, H, D, dtype=torch.float32, device=dev)
        self.rotated = w.rotated
        if self.rotated:
            # rotated basis (one per layer and KV head, shared by the sequences):
            # calibration once, then every layer's store holds the planes of (k - mu) V
            nh = w.kv_heads
            calib = torch.stack([synth.unit_calib(w, g, dev) for g in range(w.layers * nh)]).contiguous()
            self.kmean, self.kV, lam = B.fathom_calibrate_klt(calib)
            del calib
        for l in range(L):
            units = w.layer_units(l)
            keys = torch.stack([synth.unit_keys(w, u, dev) for u in units]).to(torch.bfloat16)
            if self.rotated:
                g0 = l * nh
                rk = B.fathom_rotate_keys(self.shape, keys, nh, self.kmean[g0:g0 + nh], self.kV[g0:g0 + nh])
                p, s = B.fathom_quantize_pack(self.shape, rk)
                if l == 0:
                    self.rkeys = rk                    # the rotated keys layer 0's store was coded from
                del rk
                self.var[l] = lam[g0:g0 + nh].repeat(H // nh, 1)    # unit i of the layer: head i % nh
            else:
                p, s = B.fathom_quantize_pack(self.shape, keys)
                calib = torch.stack([synth.unit_calib(w, u, dev) for u in units])
                _, self.var[l] = B.fathom_calibrate(calib)
            self.planes[l].copy_(p)
            self.scales[l].copy_(s)
            self.krows[l].copy_(keys)
            del keys, p, s
            vals = torch.stack([synth.unit_values(w, u, dev) for u in units]).to(torch.bfloat16)
            self.vrows[l].copy_(vals)
            del vals
        torch.cuda.synchronize()
        log(f"[bench] store built in {time.time() - t0:.1f}s "
            f"({'pinned host' if self.host else 'HBM'}: store {self.planes.numel() * 8 / 2**30:.2f} GiB "
            f"+ {self.scales.numel() * 2 / 2**30:.2f} GiB, rows {2 * self.krows.numel() * 2 / 2**30:.2f} GiB)")
        # queries of every step and layer (device) and their pinned host copy
        self.Q = torch.stack([torch.stack([torch.stack([synth.unit_query(w, u, dev, step=s + 1) for u in w.layer_units(l)])
                                           for l in range(L)]) for s in range(steps_total)]).contiguous()
        self.Qh = torch.empty(self.Q.shape, dtype=self.Q.dtype, pin_memory=True)
        self.Qh.copy_(self.Q)
        # per-layer budgets B_l when the workload has them (and no flat override), else flat
        self.per_layer = w.per_layer and budget <= 0
        lb = [w.budgets[l % len(w.budgets)] if self.per_layer else budget for l in range(L)]
        self.budgets = lb
        self.budget_t = torch.tensor([[b] * H for b in lb], dtype=torch.int32, device=dev)
        self.qrot = torch.empty(L, H, self.G, D, dtype=torch.float32, device=dev) if self.rotated else None
        bmax = 128 if fixed else max(lb)
        self.stage_w = max(2, min(bmax, 4 * D) * nb + (min(bmax, 4 * D) * nb) % 2)
        self.stage_s = max(8, (min(bmax, D) * nb + 7) // 8 * 8)
        self.stage_p = torch.zeros(H, self.stage_w, dtype=torch.int64, device=dev)
        self.stage_sc = torch.zeros(H, self.stage_s, dtype=torch.int16, device=dev)
        self.ws = B.alloc_workspace(self.shape, B.WS_SCAN_TOPK)
        self.aws = B.alloc_workspace(self.shape, B.WS_SPARSE_ATTN)
        self.path = path if self.host else "hbm"
        n_groups = max(1, min(groups, H))
        edges = [round(i * H / n_groups) for i in range(n_groups + 1)]
        self.groups = [(edges[i], edges[i + 1]) for i in range(n_groups) if edges[i + 1] > edges[i]]
        gsize = self.groups[0][1] - self.groups[0][0]
        assert all(b - a == gsize for a, b in self.groups), "unit groups must be equal"
        self.gshape = B.make_shape(gsize, self.n, self.D, self.G, self.k, w.n_sink, w.n_recent)
        self.gws = B.alloc_workspace(self.gshape, B.WS_SCAN_TOPK)
        self.gstream = torch.cuda.Stream()
        self.gev = [torch.cuda.Event() for _ in self.groups]
        self.depth = torch.empty(H, D, dtype=torch.uint8, device=dev)
        self.theta = torch.empty(H, dtype=torch.float64, device=dev)
        self.runs = torch.empty(H, D, 6, dtype=torch.int32, device=dev)
        self.idx = torch.empty(H, self.G, self.k, dtype=torch.int32, device=dev)
        self.sel = torch.empty(H, self.G, self.k, dtype=torch.float32, device=dev)
        self.out = torch.empty(L, H, self.G, D, dtype=torch.float32, device=dev)
        self.outh = torch.empty(L, H, self.G, D, dtype=torch.float32, pin_memory=True)
        self.qcur = torch.empty(L, H, self.G, D, dtype=torch.float32, device=dev)

    def layer(self, l, q, ev=None):
        """One layer of the decode step; ev = optional (start, end) events around the
        dominant stage (host regime: the gather, or the fused scan; HBM regime: the scan).
        A rotated store is planned and scanned with the rotated queries q V; the exact
        attention takes the original q."""
        B = self.B
        qa = q
        if self.rotated:
            nh = self.w.kv_heads
            q = B.fathom_rotate_query(self.shape, qa, nh, self.kV[l * nh:(l + 1) * nh], out=self.qrot[l])
        if self.fixed:
            B.fathom_plan_fixed(self.shape, q, self.var[l], 32, 4, depth=self.depth, runs=self.runs)
        else:
            B.fathom_plan(self.shape, q, self.var[l], self.budget_t[l], depth=self.depth, theta=self.theta,
                          runs=self.runs, want_theta=self.want_theta)
        if self.host and self.path == "pipelined":
            self._gather_scan_pipelined(l, q, ev)
        elif self.host and self.path == "staged":
            if ev:
                ev[0].record()
            B.fathom_gather(self.shape, self.planes[l], self.scales[l], self.runs, self.stage_p, self.stage_sc)
            if ev:
                ev[1].record()
            B.fathom_scan_topk(self.shape, self.stage_p, self.stage_sc, self.runs, q, self.ws,
                               source=B.SRC_STAGING, topk_idx=self.idx, topk_score=self.sel)
        else:
            # HBM regime, or the fused host path: the scan stages the planned runs
            # straight from the store (pinned host memory) into shared memory
            if ev:
                ev[0].record()
            B.fathom_scan_topk(self.shape, self.planes[l], self.scales[l], self.runs, q, self.ws,
                               topk_idx=self.idx, topk_score=self.sel)
            if ev:
                ev[1].record()
        B.fathom_sparse_attn(self.shape, self.krows[l], self.vrows[l], qa, self.idx, self.aws, out=self.out[l])

    def _gather_scan_pipelined(self, l, q, ev=None):
        """Gathers of unit groups on a second stream, each group's scan on the main stream
        as soon as its runs have landed in HBM staging: the link stays busy while the SMs scan."""
        B = self.B
        main = torch.cuda.current_stream()
        gs = self.gstream
        plan_done = torch.cuda.Event()
        plan_done.record(main)             # also orders this layer's gathers after the last layer's scans
        gs.wait_event(plan_done)
        n_g = len(self.groups)
        if ev:
            ev[0].record(gs)
        for g, (a, b) in enumerate(self.groups):
            with torch.cuda.stream(gs):
                B.fathom_gather(self.gshape, self.planes[l, a:b], self.scales[l, a:b], self.runs[a:b],
                                self.stage_p[a:b], self.stage_sc[a:b])
                if ev and g == n_g - 1:
                    ev[1].record(gs)
                self.gev[g].record(gs)
            main.wait_event(self.gev[g])
            B.fathom_scan_topk(self.gshape, self.stage_p[a:b], self.stage_sc[a:b], self.runs[a:b], q[a:b],
                               self.gws, source=B.SRC_STAGING, topk_idx=self.idx[a:b], topk_score=self.sel[a:b])

    def layer_stages(self, l, q):
        """One layer with CUDA events between the calls: per-stage milliseconds (the
        pipelined path reports its overlapped gather + scan as one stage)."""
        B = self.B
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        qa = q
        ev[0].record()
        if self.rotated:
            nh = self.w.kv_heads
            q = B.fathom_rotate_query(self.shape, qa, nh, self.kV[l * nh:(l + 1) * nh], out=self.qrot[l])
        if self.fixed:
            B.fathom_plan_fixed(self.shape, q, self.var[l], 32, 4, depth=self.depth, runs=self.runs)
        else:
            B.fathom_plan(self.shape, q, self.var[l], self.budget_t[l], depth=self.depth, theta=self.theta,
                          runs=self.runs, want_theta=self.want_theta)
        ev[1].record()
        if self.host and self.path == "staged":
            B.fathom_gather(self.shape, self.planes[l], self.scales[l], self.runs, self.stage_p, self.stage_sc)
            ev[2].record()
            B.fathom_scan_topk(self.shape, self.stage_p, self.stage_sc, self.runs, q, self.ws,
                               source=B.SRC_STAGING, topk_idx=self.idx, topk_score=self.sel)
        elif self.host and self.path == "pipelined":
            ev[2].record()
            self._gather_scan_pipelined(l, q)
        else:
            ev[2].record()
            B.fathom_scan_topk(self.shape, self.planes[l], self.scales[l], self.runs, q, self.ws,
                               topk_idx=self.idx, topk_score=self.sel)
        ev[3].record()
        B.fathom_sparse_attn(self.shape, self.krows[l], self.vrows[l], qa, self.idx, self.aws, out=self.out[l])
        ev[4].record()
        return ev

    def capture(self, evs):
        """One decode step (all layers) as a CUDA graph reading the queries from
        self.qcur; evs[l] = events (recorded inside the graph) around layer l's
        dominant stage."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):          # warm the calls on the capture stream's side
            for l in range(self.L):
                self.layer(l, self.qcur[l])
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for l in range(self.L):
                self.layer(l, self.qcur[l], evs[l] if evs else None)
        torch.cuda.synchronize()
        return g

    def step(self, s, evs=None):
        for l in range(self.L):
            self.layer(l, self.Q[s, l], evs[l] if evs else None)

    def step_e2e(self, s):
        """The same step through the public calls with host buffers: the step's
        queries come from pinned host memory and the attention outputs go back."""
        self.qcur.copy_(self.Qh[s], non_blocking=True)
        for l in range(self.L):
            self.layer(l, self.qcur[l])
        self.outh.copy_(self.out, non_blocking=True)

    def planned_bytes(self):
        """Scanned bytes of the current plan per layer (code planes + active scales), summed over units."""
        d = self.depth.to(torch.int64)
        return int(d.sum().item()) * self.nb * 8 + int((d > 0).sum().item()) * self.nb * 2


def measure_link_peak():
    """Pinned host -> device copy bandwidth (copy engine), best of 10 over 1 GiB."""
    sz = 1 << 30
    h = torch.empty(sz, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(sz, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    best = 1e9
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / 1e3)
    del h, d
    return sz / best / 1e9


def measure_sm_read_peak(st):
    """Host-link read rate of SM loads (not the copy engine): fathom_gather of a plan with
    every channel at depth 4 copies layer 0's whole pinned store (68 B per token and unit)
    into HBM with 16-byte loads from every SM; best of 5."""
    B = st.B
    H, D, nb = st.H, st.D, st.nb
    q = st.Q[0, 0]
    depth, runs = B.fathom_plan_fixed(st.shape, q, st.var[0], D, 4)
    sp = torch.empty(H, 4 * D * nb, dtype=torch.int64, device="cuda")
    ss = torch.empty(H, D * nb + (-(D * nb)) % 8, dtype=torch.int16, device="cuda")
    nbytes = H * (4 * D * nb * 8 + D * nb * 2)
    for _ in range(2):
        B.fathom_gather(st.shape, st.planes[0], st.scales[0], runs, sp, ss)
    torch.cuda.synchronize()
    best = 1e9
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        B.fathom_gather(st.shape, st.planes[0], st.scales[0], runs, sp, ss)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / 1e3)
    del sp, ss
    return nbytes / best / 1e9


# Thread instructions the first-pass scan kernel issues per scored token, from the
# ncu capture of one HBM-resident host_1m layer (8 units x 2^20 tokens, B = 48) of
# the current kernel; the bench multiplies it by the tokens a call scores to
# estimate how close the HBM-resident scan runs to the instruction-issue bound.
SCAN_PROFILE = {"thread_instructions_per_token": 71.59e6 * 32 / (8 << 20),
                "dram_bytes_per_layer": 56.98e6 + 0.87e6,
                "source": "profiles/scan_kernel_host1m_hbm.md"}


def measure_hbm_scan(st, args, peaks, sm_mhz):
    """The scan + top-k call on layer 0's store copied into HBM (the HBM-resident
    regime), with each timed step's plan; L2 (129 MB) is flushed by a 256 MiB write
    before every call, and CUDA events bracket the call on its stream."""
    B = st.B
    planes = st.planes[0].to("cuda")
    scales = st.scales[0].to("cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    times, nbytes = [], []
    for i in range(args.warmup + args.steps):
        q = st.Q[i, 0]
        if st.fixed:
            B.fathom_plan_fixed(st.shape, q, st.var[0], 32, 4, depth=st.depth, runs=st.runs)
        else:
            B.fathom_plan(st.shape, q, st.var[0], st.budget_t[0], depth=st.depth, runs=st.runs, want_theta=False)
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        B.fathom_scan_topk(st.shape, planes, scales, st.runs, q, st.ws, topk_idx=st.idx, topk_score=st.sel)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
            nbytes.append(st.planned_bytes())
    del planes, scales, flush
    t = statistics.mean(times)
    gbs = statistics.mean(nbytes) / t / 1e9
    hbm = peaks["hbm_gbs"]
    res = {"us": t * 1e6, "gbs": gbs, "peak_gbs": hbm, "frac": gbs / hbm,
           "scanned_bytes": statistics.mean(nbytes), "calls": len(times),
           "traffic": SCAN_PROFILE["dram_bytes_per_layer"],
           "note": "fathom_scan_topk (first-pass scan, merge, exact second pass, second merge) on layer 0's "
                   "store copied to HBM, the plan of each timed step's queries, L2 flushed before each call; "
                   "traffic = DRAM read + write bytes of the first-pass scan kernel on this layer "
                   f"({SCAN_PROFILE['source']})"}
    ipt = SCAN_PROFILE["thread_instructions_per_token"]
    if ipt:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        mhz = sm_mhz or 2070.0
        tokens = st.H * st.n
        res["issue_bound_frac"] = ipt * tokens / 32.0 / (sms * 4 * mhz * 1e6 * t)
        res["issue_note"] = (f"{ipt:.0f} thread instructions per token (profiled) x {tokens} tokens / 32 = warp "
                             f"instructions, over {sms} SMs x 4 issue slots x {mhz:.0f} MHz x the call's time")
    return res


def measure_fixed_plan(st, args):
    """The byte-equivalent 136-bit comparison (32 channels at depth 4, the same kernels),
    timed as the main step: one graph replay per step, each with its own queries."""
    st.fixed = True
    try:
        graph = st.capture(None)
        gw = max(args.warmup, 10)
        for i in range(gw):
            st.qcur.copy_(st.Q[i], non_blocking=True)
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(args.steps):
            st.qcur.copy_(st.Q[gw + i], non_blocking=True)
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        us_layer = e0.elapsed_time(e1) * 1e3 / (args.steps * st.L)
        st.layer(0, st.Q[0, 0])
        torch.cuda.synchronize()
        nbytes = st.planned_bytes()
        del graph
    finally:
        st.fixed = False
    return {"us_per_layer": us_layer, "scanned_bytes_per_layer": nbytes}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return json.load(open(p)), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ---------------------------------------------------------------- CPU oracle baseline
def unit_budget(w: synth.Workload, budget: int, unit: int) -> int:
    """The unit's code-bit budget: the flat budget, or its layer's B_l (budget <= 0)."""
    if w.per_layer and budget <= 0:
        return w.budgets[((unit // w.kv_heads) % w.layers) % len(w.budgets)]
    return budget


def _oracle_inputs(w: synth.Workload, budget: int, unit: int) -> dict:
    """One unit's inputs to the oracle's decode step, with its store built (the
    store build is not part of the step and is not timed)."""
    from oracle import oracle as O
    O.build()
    keys = synth.unit_keys(w, unit, "cpu").to(torch.bfloat16)
    k32 = keys.float().numpy()
    kb = keys.view(torch.int16).numpy().view(np.uint16)
    vb = synth.unit_values(w, unit, "cpu").to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q = synth.unit_query(w, unit, "cpu", step=1).numpy()
    calib = synth.unit_calib(w, unit, "cpu").numpy()
    V = None
    if w.rotated:
        mean, _, cov = O.calibrate(calib, with_cov=True)
        lam, V = O.eigh(cov)
        var = lam.astype(np.float32)
        k32 = O.rotate(k32, mean, V)
    else:
        _, var = O.calibrate(calib)
        var = var.astype(np.float32)
    P, S, _ = O.quantize_pack(k32)
    return {"kb": kb, "vb": vb, "q": q, "V": V, "var": var, "P": P, "S": S,
            "budget": unit_budget(w, budget, unit)}


def _oracle_step(w: synth.Workload, inp: dict) -> float:
    """The oracle's whole per-unit decode step (query rotation for a rotated
    store, plan, gather, scores, selection, attention); returns seconds."""
    from oracle import oracle as O
    n = w.n
    t0 = time.perf_counter()
    qs = O.rotate_query(inp["q"], inp["V"]).astype(np.float32) if w.rotated else inp["q"]
    depth, theta, _ = O.plan(qs, inp["var"], inp["budget"])
    runs = O.runs(depth, n)
    if w.regime == "host":
        nb = (n + 63) // 64
        sp, ss = O.gather(runs, inp["P"], inp["S"], int(depth.sum()) * nb, int((depth > 0).sum()) * nb)
        s = O.scores_staged(runs, sp, ss, depth, qs, n)
    else:
        s = O.scores(inp["P"][None], inp["S"][None], depth[None], qs[None], n)[0]
    idx, _ = O.select(s, w.k, w.n_sink, w.n_recent)
    O.attention(inp["kb"], inp["vb"], inp["q"], idx)
    return time.perf_counter() - t0


def oracle_layer_sample(w: synth.Workload, budget: int, unit: int):
    """Time the CPU oracle on one unit of the workload; returns seconds."""
    return _oracle_step(w, _oracle_inputs(w, budget, unit))


def cpu_baseline(w, budget, reps=1):
    secs = [oracle_layer_sample(w, budget, u) for u in w.layer_units(0)[:reps]]
    per_unit = statistics.mean(secs)
    us_layer = per_unit * w.units_per_layer() * 1e6
    return {"value": us_layer, "unit": "µs/layer", "cores": 1, "kind": "oracle",
            "sample": f"{reps} unit(s) of layer 0 at n={w.n} (plan, gather, scores, top-k, attention; "
                      f"single-threaded C), scaled x{w.units_per_layer()} units per layer"}


def _parallel_worker(w: synth.Workload, budget: int, unit: int, barrier, wait_s: float, results):
    """One worker process of the all-cores baseline: build the unit's inputs,
    wait for the other workers, then time the unit's step (monotonic clock,
    comparable across the processes of one host).  Puts (unit, t0, t1) or
    (unit, error) on `results`."""
    try:
        torch.set_num_threads(1)
        inp = _oracle_inputs(w, budget, unit)
        barrier.wait(timeout=wait_s)
        t0 = time.monotonic()
        _oracle_step(w, inp)
        results.put((unit, t0, time.monotonic()))
    except BaseException as exc:   # the parent reports it; never hang the barrier's other parties
        try:
            barrier.abort()
        finally:
            results.put((unit, repr(exc)[:200]))


def host_cores() -> int:
    """Cores this process may run on (its affinity set)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline_parallel(w: synth.Workload, budget: int, max_workers: int = 0, mem_bytes: int = 8 << 30,
                          wait_s: float = 600.0) -> dict:
    """The oracle on several units of layer 0 at once, one single-threaded process per
    unit ("spawn" processes: this process already holds a CUDA context).  Workers are
    limited by the host's cores, the layer's units and a host-memory budget for their
    inputs (about 14 bytes per token and channel).  The layer's time is the wall time
    of one round (first start to last end, after a barrier) times the rounds a layer
    needs on that many workers.  A worker that fails or does not report within
    2 * wait_s is terminated and the call raises."""
    import math
    import multiprocessing as mp
    import queue as queue_mod
    per_unit = 14 * w.n * w.D
    P = min(host_cores(), w.units_per_layer(), max(1, mem_bytes // per_unit))
    if max_workers:
        P = min(P, max_workers)
    P = max(1, P)
    units = w.layer_units(0)[:P]
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(P), ctx.Queue()
    procs = [ctx.Process(target=_parallel_worker, args=(w, budget, u, barrier, wait_s, results), daemon=True)
             for u in units]
    spans, errors = [], []
    try:
        for pr in procs:
            pr.start()
        deadline = time.monotonic() + 2 * wait_s
        while len(spans) + len(errors) < P:
            try:
                r = results.get(timeout=2.0)
            except queue_mod.Empty:
                dead = [pr.exitcode for pr in procs if not pr.is_alive() and pr.exitcode not in (0, None)]
                if dead:
                    raise RuntimeError(f"all-cores baseline: a worker exited with code {dead[0]}")
                if time.monotonic() > deadline:
                    raise TimeoutError(f"all-cores baseline: {P - len(spans) - len(errors)} worker(s) "
                                       "did not report")
                continue
            (spans if len(r) == 3 else errors).append(r)
    finally:
        for pr in procs:
            pr.join(timeout=10)
            if pr.is_alive():
                pr.terminate()
                pr.join(timeout=10)
    if errors:
        raise RuntimeError(f"all-cores baseline: worker error {errors[0]}")
    wall = max(t1 for _, _, t1 in spans) - min(t0 for _, t0, _ in spans)
    rounds = math.ceil(w.units_per_layer() / P)
    return {"value": wall * rounds * 1e6, "unit": "µs/layer", "cores": P, "kind": "oracle",
            "sample": f"{P} unit(s) of layer 0 at n={w.n} in {P} single-threaded processes at once "
                      f"(wall time of the round), x{rounds} rounds for the layer's "
                      f"{w.units_per_layer()} units; {host_cores()} cores available"}


# ---------------------------------------------------------------- main
def workload_config(w: synth.Workload, args) -> dict:
    """The JSON line's config (the same for both arms)."""
    per_layer = w.per_layer and args.budget <= 0
    budgets = [w.budgets[l % len(w.budgets)] if per_layer else args.budget for l in range(w.layers)]
    path = args.path if w.regime == "host" else "hbm"
    return {"workload": w.name, "n": w.n, "layers": w.layers, "kv_heads": w.kv_heads, "sessions_per_gpu": w.seqs,
            "G": w.G, "D": w.D, "k": w.k, "n_sink": w.n_sink, "n_recent": w.n_recent,
            "budget": ("fixed 32ch x 4 planes" if args.fixed else
                       f"per layer {budgets}" if per_layer else args.budget),
            "basis": "rotated (KLT per layer and KV head)" if w.rotated else "channels",
            "regime": w.regime, "path": path,
            "unit_groups": args.groups if path == "pipelined" else 1,
            "l2": l2_note(w)}


L2_BYTES = 129 << 20      # GB300 L2
# Graph replays before the timed region.  On a host-resident store the first
# replays run slower (up to 1.4x over the first ten or so, in every run) while
# the pinned pages' translations warm up; a decode loop runs in the steady state
# that follows.
GRAPH_WARMUP = 40


def l2_note(w: synth.Workload) -> str:
    """Whether the step's inputs exceed L2 (the timing rule: inputs larger than L2,
    or an L2 flush between timed steps; this bench never flushes)."""
    store = w.units * w.n * (w.D // 2 + w.D // 32)      # 4 plane bits + a 16-bit scale per 64 tokens
    rows = w.units * w.n * w.D * 2 * 2                   # bf16 K and V rows
    mb = (store + rows) / 2**20
    if store + rows > L2_BYTES:
        return f"inputs larger than L2 (store and rows of all layers: {mb:.0f} MiB > 129 MiB)"
    return f"inputs fit in L2 ({mb:.1f} MiB): L2-resident, latency-bound; no HBM roofline claim"


def run_reference(args, w, rank, world):
    """The CPU oracle on the same workload, as the reference arm.  One step is one
    (layer, KV head) unit's decode step, which is what is timed: ms_per_step is that
    unit's time, and value scales it to a layer (x units per layer) so that it
    reads in the same unit as the GPU arm's value."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_layer_sample(w, args.budget, w.layer_units(0)[0])
    secs = []
    units = w.layer_units(0)
    for s in range(args.steps):
        secs.append(oracle_layer_sample(w, args.budget, units[s % len(units)]))
    per_unit = statistics.mean(secs)
    us_layer = per_unit * w.units_per_layer() * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": us_layer, "unit": "µs/layer",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_unit * 1e3,
            "step": f"one unit (one KV head of one layer) at n={w.n}; value = the unit's time x "
                    f"{w.units_per_layer()} units per layer",
            "unit_step_ms_min_median_max": [min(secs) * 1e3, statistics.median(secs) * 1e3, max(secs) * 1e3],
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Qwen3-8B-shaped keys/queries/values)",
            "config": workload_config(w, args),
            "cpu_baseline": {"value": us_layer, "unit": "µs/layer", "cores": 1, "kind": "oracle",
                             "sample": f"one unit per step at n={w.n}, scaled x{w.units_per_layer()} units per layer"},
            "e2e": {"value": us_layer, "unit": "µs/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def spawn_ranks(n):
    """`--gpus N` without a launcher: start N copies of this command as ranks
    0..N-1 of one job on this node (RANK, LOCAL_RANK, WORLD_SIZE and a free
    MASTER_PORT on 127.0.0.1 in their environment), pass rank 0's output
    through, and return the largest exit code."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    procs = []
    for r in range(n):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        out = None if r == 0 else subprocess.DEVNULL
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__), *sys.argv[1:]], env=env,
                                      stdout=out))
    rcs = [p.wait() for p in procs]
    return max(abs(rc) for rc in rcs)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="host_1m", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--budget", type=int, default=None,
                    help="flat code-bit budget (default: 48, or the per-layer budgets of a workload that has them)")
    ap.add_argument("--fixed", action="store_true", help="the 136-bit fixed-depth comparison plan")
    ap.add_argument("--path", default="fused", choices=["fused", "staged", "pipelined"],
                    help="host regime: the scan reads the pinned store directly (default), gather then "
                         "scan, or gathers overlapped with scans")
    ap.add_argument("--groups", type=int, default=4, help="unit groups of the pipelined path")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of a CUDA graph per step")
    ap.add_argument("--impl", default="fathom", choices=["fathom", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (0: workload's)")
    ap.add_argument("--regime", default="", choices=["", "hbm", "host"],
                    help="override where the store and rows live (default: the workload's)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fidelity", action="store_true", help="skip the (untimed) fidelity measurement")
    ap.add_argument("--plan-theta", action="store_true",
                    help="have the plan also write theta (the decode step needs only the depths and runs)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the HBM-resident scan and 136-bit comparison measurements")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_ranks(args.gpus))
    if int(os.environ.get("WORLD_SIZE", "1")) != args.gpus:
        log(f"[bench] --gpus {args.gpus} but WORLD_SIZE={os.environ.get('WORLD_SIZE')}: launch one rank per GPU")
        sys.exit(2)
    rank, world = dist_setup(args.gpus)
    w = synth.WORKLOADS[args.workload]
    if args.budget is None:
        args.budget = 0 if w.per_layer else 48
    if args.layers:
        w = synth.shrink(w, layers=args.layers)
    if args.regime:
        w = synth.shrink(w, regime=args.regime)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    from bit_plane_kv_gb300 import binding as B
    import __graft_entry__
    __graft_entry__.build()
    # queries: warm-up, timed, e2e, graph warm-up and 50 spread steps, all distinct
    total_steps = args.warmup + 2 * args.steps + max(args.warmup, GRAPH_WARMUP) + 50
    st = Setup(w, args.budget, rank, total_steps, args.fixed, args.path, args.groups, args.plan_theta)
    link_gbs = measure_link_peak() if st.host else None
    sm_link_gbs = measure_sm_read_peak(st) if st.host else None
    link_src = "measured in this run: pinned host->device copy, 1 GiB, best of 10"
    if st.host and sm_link_gbs > link_gbs:
        link_gbs, link_src = sm_link_gbs, "measured in this run: SM loads of the whole pinned store (fathom_gather), best of 5"
    peaks, peak_src = measured_peaks()

    # warm-up
    for s in range(args.warmup):
        st.step(s)
    torch.cuda.synchronize()
    plan_bytes = [0] * st.L
    active = [0.0] * st.L                 # mean active channels (t_j > 0) per unit, per layer
    for l in range(st.L):
        st.layer(l, st.Q[0, l])
        torch.cuda.synchronize()
        plan_bytes[l] = st.planned_bytes()
        active[l] = float((st.depth > 0).sum().item()) / st.H

    # CPU time to issue one eager step (the Python binding's per-call cost)
    torch.cuda.synchronize()
    c0 = time.perf_counter()
    st.step(0)
    issue_s = time.perf_counter() - c0
    torch.cuda.synchronize()

    # timed region: K steps, each one replay of the step's CUDA graph (queries
    # copied into the graph's input buffer first), with events captured around
    # the dominant stage of every layer
    use_graph = not args.eager
    try:
        gevs = [(torch.cuda.Event(enable_timing=True, external=True),
                 torch.cuda.Event(enable_timing=True, external=True)) for _ in range(st.L)] if use_graph else None
        graph = st.capture(gevs) if use_graph else None
    except Exception as exc:               # no graph capture: time the eager step
        log(f"[bench] CUDA graph capture unavailable ({exc}); timing eager launches")
        use_graph, graph = False, None
    clocks = ClockSampler()
    clocks.start()                              # running (first sample taken) before the timed region
    # graph warm-up: the first replays upload the graph, and a host-resident store needs
    # several steps with different queries (different planned channels) before its reads
    # reach their steady rate, as in a decode loop: at least GRAPH_WARMUP replays, each with its own
    # queries (none of them used by the timed steps)
    graph_warmup = max(args.warmup, GRAPH_WARMUP) if use_graph else 0
    q_gw = args.warmup + 2 * args.steps         # first query index reserved for the graph warm-up
    if use_graph:
        for s in range(graph_warmup):
            st.qcur.copy_(st.Q[q_gw + s], non_blocking=True)
            graph.replay()
        torch.cuda.synchronize()
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(st.L)]
           for _ in range(args.steps)]
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kern = []
    t_start.record()
    step_ev[0].record()
    for s in range(args.steps):
        if use_graph:
            st.qcur.copy_(st.Q[args.warmup + s], non_blocking=True)
            graph.replay()
        else:
            st.step(args.warmup + s, evs[s])
        step_ev[s + 1].record()
    t_end.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    clk = clocks.stop(torch.cuda.current_device(), window=(wall0, wall1))
    elapsed = t_start.elapsed_time(t_end) / 1e3
    step_ms = [step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps)]
    log("[bench] step ms: " + " ".join(f"{x:.3f}" for x in step_ms))
    elapsed = max_over_ranks(elapsed, world)
    if use_graph:
        # the captured events hold the last replay's stage times; one more replay per step for the average
        for s in range(args.steps):
            st.qcur.copy_(st.Q[args.warmup + s], non_blocking=True)
            graph.replay()
            torch.cuda.synchronize()
            kern += [a.elapsed_time(b) / 1e3 for a, b in gevs]
    else:
        kern = [e[0].elapsed_time(e[1]) / 1e3 for row in evs for e in row]
    kern_avg = statistics.mean(kern)

    # end to end through the public calls with host buffers, on the host clock: each
    # step issues its query copy, every layer's calls and the output copy, and waits
    # for the output (a decode loop reads it before the next step)
    barrier(world)
    torch.cuda.synchronize()
    e2e_steps = []
    for s in range(args.steps):
        h0 = time.perf_counter()
        st.step_e2e(args.warmup + args.steps + s)
        torch.cuda.current_stream().synchronize()
        e2e_steps.append(time.perf_counter() - h0)
    e2e_elapsed = max_over_ranks(sum(e2e_steps), world)

    # per-step spread over more steps than the timed region (graph replays, each with
    # its own queries; events between replays), reported beside the timed value
    spread_ms = []
    if use_graph:
        n_spread = 50
        sp_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_spread + 1)]
        q_sp = args.warmup + 2 * args.steps + graph_warmup
        sp_ev[0].record()
        for i in range(n_spread):
            st.qcur.copy_(st.Q[q_sp + i], non_blocking=True)
            graph.replay()
            sp_ev[i + 1].record()
        torch.cuda.synchronize()
        spread_ms = sorted(sp_ev[i].elapsed_time(sp_ev[i + 1]) for i in range(n_spread))

    # decode-time append: coding the block of a new token into the store (the step before
    # the scan in a decode loop); timed on layer 0's store for its last block, which codes
    # the same values again, as a graph of `steps` appends
    append_us = None
    try:
        B = st.B
        blk, cnt = (st.n - 1) // 64, (st.n - 1) % 64 + 1
        keys_l0 = st.rkeys if st.rotated else st.krows[0]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            B.fathom_append_block(st.shape, keys_l0, blk, cnt, st.planes[0], st.scales[0])
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        ag = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ag):
            for _ in range(args.steps):
                B.fathom_append_block(st.shape, keys_l0, blk, cnt, st.planes[0], st.scales[0])
        ag.replay()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        ag.replay()
        a1.record()
        torch.cuda.synchronize()
        append_us = a0.elapsed_time(a1) * 1e3 / args.steps
    except Exception as exc:   # reported as missing, never as a number
        log(f"[bench] append timing unavailable: {exc}")

    # the HBM-resident scan and the 136-bit comparison (host-resident runs)
    hbm_scan, fixed136 = None, None
    if st.host and not args.no_extras:
        try:
            hbm_scan = measure_hbm_scan(st, args, peaks, clk.get("sm_mhz"))
            log(f"[bench] HBM-resident scan: {hbm_scan}")
        except Exception as exc:   # reported as missing, never as a number
            log(f"[bench] HBM-resident scan unavailable: {exc}")
            hbm_scan = {"error": str(exc)[:200]}
        if not st.fixed and st.path == "fused":
            try:
                fixed136 = measure_fixed_plan(st, args)
                log(f"[bench] 136-bit plan: {fixed136}")
            except Exception as exc:   # reported as missing, never as a number
                log(f"[bench] 136-bit plan unavailable: {exc}")
                fixed136 = {"error": str(exc)[:200]}

    # per-stage breakdown (separate pass, events between the calls)
    stage_ev = []
    for s in range(args.steps):
        for l in range(st.L):
            stage_ev.append(st.layer_stages(l, st.Q[args.warmup + s, l]))
    torch.cuda.synchronize()
    names = ["plan", "gather", "scan_topk", "sparse_attn"]
    stages = {nm: statistics.mean(e[i].elapsed_time(e[i + 1]) * 1e3 for e in stage_ev) for i, nm in enumerate(names)}
    log("[bench] per-layer stages (µs): " + ", ".join(f"{k} {v:.1f}" for k, v in stages.items()))

    # rotated workloads: the calibration-free basis from the sessions' own keys
    # (one layer of the workload, and one layer of 8 KV heads at 100k tokens)
    klt_online = None
    if st.rotated:
        try:
            B = st.B

            def time_online(shape, rows, reps=3):
                ws = B.alloc_workspace(shape, B.WS_KLT_ONLINE)
                m = torch.empty(shape.units, shape.D, dtype=torch.float64, device="cuda")
                V = torch.empty(shape.units, shape.D, shape.D, dtype=torch.float64, device="cuda")
                lam = torch.empty(shape.units, shape.D, dtype=torch.float32, device="cuda")
                for _ in range(2):
                    B.fathom_klt_online(shape, rows, ws, m, V, lam)
                torch.cuda.synchronize()
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record()
                for _ in range(reps):
                    B.fathom_klt_online(shape, rows, ws, m, V, lam)
                a1.record()
                torch.cuda.synchronize()
                return a0.elapsed_time(a1) * 1e3 / reps

            us_layer = time_online(st.shape, st.krows[0])
            units8 = st.w.layer_units(0)[:8]
            rows100k = torch.stack([synth.unit_keys(st.w, u, "cuda", n=100000) for u in units8]).to(torch.bfloat16)
            us_100k = time_online(B.make_shape(8, 100000, st.D, st.G, 1, 0, 0), rows100k)
            del rows100k
            klt_online = {"us_per_layer": us_layer, "layer_units": st.H, "layer_tokens": st.n,
                          "us_8_heads_100k_tokens": us_100k,
                          "note": "fathom_klt_online (mean, covariance, fp32 Jacobi) on each unit's own keys, "
                                  "CUDA events, mean of 3 calls after 2 warm-up calls"}
            log(f"[bench] online basis: {klt_online}")
        except Exception as exc:   # reported as missing, never as a number
            log(f"[bench] online basis timing unavailable: {exc}")
            klt_online = {"error": str(exc)[:200]}

    # fidelity of the timed path (untimed): layer 0 at the last timed step's query,
    # against dense attention and against attention over the exact top-k
    fidelity = None
    if not args.no_fidelity:
        try:
            from bit_plane_kv_gb300 import fidelity as FID
            q0 = st.Q[args.warmup + args.steps - 1, 0].contiguous()
            st.layer(0, q0)
            res = FID.compare(st.shape, st.krows[0], st.vrows[0], q0, st.idx, st.out[0],
                              workspaces={"scan": st.ws, "attn": st.aws})
            # the same kept sets attended with keys rebuilt from the store's four planes
            # (no bf16 K rows), timed over 3 calls
            B = st.B
            qk = st.qrot[0] if st.rotated else q0
            pl_out = torch.empty_like(st.out[0])
            B.fathom_sparse_attn_planes(st.shape, st.planes[0], st.scales[0], st.vrows[0], qk, st.idx, st.aws, out=pl_out)
            torch.cuda.synchronize()
            p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            p0.record()
            for _ in range(3):
                B.fathom_sparse_attn_planes(st.shape, st.planes[0], st.scales[0], st.vrows[0], qk, st.idx, st.aws,
                                            out=pl_out)
            p1.record()
            torch.cuda.synchronize()
            dense0 = B.fathom_dense_attn(st.shape, st.krows[0], st.vrows[0], q0,
                                         B.alloc_workspace(st.shape, B.WS_DENSE_ATTN))
            rel_pl = B.fathom_rel_err(pl_out, dense0).cpu().numpy()
            rel_pl_rows = B.fathom_rel_err(pl_out, st.out[0]).cpu().numpy()
            fidelity = {
                "layer": 0, "budget": st.budgets[0] if not st.fixed else "fixed 136-bit",
                "planes_k_rel_l2_vs_dense_mean": float(rel_pl.mean()),
                "planes_k_rel_l2_vs_bf16_k_mean": float(rel_pl_rows.mean()),
                "planes_k_attn_us_per_layer": p0.elapsed_time(p1) * 1e3 / 3,
                "rel_l2_vs_dense_mean": float(res["rel_dense"].mean()),
                "rel_l2_vs_dense_max": float(res["rel_dense"].max()),
                "rel_l2_vs_exact_topk_mean": float(res["rel_exact"].mean()),
                "exact_topk_rel_l2_vs_dense_mean": float(res["exact_vs_dense"].mean()),
                "exact_topk_overlap_mean": float(res["overlap"].mean()),
                "note": "relative L2 error of the attention output per (unit, head), averaged; overlap = "
                        "fraction of the exact top-k (q . k over the bf16 rows) the scan kept; planes_k: the "
                        "kept sets attended with keys rebuilt from the store's four planes instead of bf16 K rows",
            }
            log(f"[bench] fidelity: {fidelity}")
        except Exception as exc:   # reported as missing, never as a number
            log(f"[bench] fidelity unavailable: {exc}")
            fidelity = {"error": str(exc)[:200]}

    L, H = st.L, st.H
    layer_steps = args.steps * L * world
    us_layer = elapsed * 1e6 / layer_steps         # whole job: all ranks' layer-steps
    e2e_us_layer = e2e_elapsed * 1e6 / layer_steps
    scanned = statistics.mean(plan_bytes)          # bytes scanned per layer (all units of the layer)
    bits_per_token = scanned * 8 / (H * st.n)
    scan_gbs = scanned / (elapsed / (args.steps * L)) / 1e9
    # our kernel launches per layer: plan, attention, and scan_topk's four (scan,
    # merge, exact second-pass scan, second merge), plus one gather per group
    if st.host and st.path == "pipelined":
        launches_per_layer = 2 + 5 * len(st.groups)
    elif st.host and st.path == "staged":
        launches_per_layer = 7
    else:
        launches_per_layer = 6
    launches_per_layer += 1 if st.rotated else 0     # the query rotation
    if st.host:
        link = link_gbs
        achieved = scanned / kern_avg / 1e9
        what = {"staged": ("gather_kernel", "gather launch"),
                "pipelined": ("gather_kernel", "layer's gather launches (one per unit group, back to back on "
                                               "their own stream, overlapped with the scans)"),
                "fused": ("scan_kernel", "fused scan_topk call (its scan kernel loads the runs from pinned "
                                         "host memory)")}[st.path]
        roof = {"bound": "link", "achieved": achieved, "peak": link, "unit": "GB/s", "frac": achieved / link,
                "traffic": None, "kernel": what[0],
                "traffic_note": "the runs cross the host link, not HBM: no DRAM counter measures them",
                "peak_source": link_src + " (the larger of the copy-engine and SM-load rates)",
                "note": f"host-link bytes (planned plane runs + active-channel scales) per {what[1]} / its time"}
    else:
        hbm = peaks["hbm_gbs"]
        achieved = scanned / kern_avg / 1e9
        same_as_profile = w.name == "host_1m" and args.budget == 48 and not args.fixed
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": SCAN_PROFILE["dram_bytes_per_layer"] if same_as_profile else None,
                "kernel": "scan_kernel",
                "traffic_note": (f"DRAM read + write bytes of the first-pass scan kernel on one layer of this "
                                 f"workload ({SCAN_PROFILE['source']})" if same_as_profile else
                                 "no ncu capture of this workload's scan layer"),
                "peak_source": f"{peak_src} HBM copy peak (MEASURED_PEAKS.json hbm_gbs)",
                "binding_resource": f"instruction issue ({SCAN_PROFILE['source']})",
                "note": "scanned bytes per layer / the scan_topk call's time (scan + merge kernels); the HBM "
                        "roofline is the denominator the target is stated against, not the scan's bound"}
    line = {
        "metric": METRIC, "value": us_layer, "unit": "µs/layer", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp32 (u64 bit planes, fp16 scales, bf16 rows)",
        "data": "synthetic (seeded Qwen3-8B-shaped keys/queries/values, no trained weights)",
        "config": workload_config(w, args),
        "scan_gbs": scan_gbs,
        "scanned_bytes_per_layer": scanned,
        "scanned_bits_per_token": bits_per_token,
        "active_channels_per_unit": statistics.mean(active),
        "roofline": roof,
        "e2e": {"value": e2e_us_layer, "unit": "µs/layer",
                "h2d_bytes_per_step": int(st.Q[0].numel() * 4), "d2h_bytes_per_step": int(st.out.numel() * 4),
                "how": "host wall clock (perf_counter) per step around the query copy from pinned host memory, "
                       "every layer's C-ABI calls (eager, through the Python binding) and the output copy back, "
                       "ending at the stream's synchronisation"},
        "gpu_launches": launches_per_layer * L * args.steps,
        "stages_us_per_layer": stages,
        "append_us_per_layer": append_us,
        "fidelity": fidelity,
        "klt_online": klt_online,
        "timing": "one CUDA graph replay per step" if use_graph else "eager launches",
        "graph_warmup_replays": graph_warmup,
        "step_ms_min_median_max": [min(step_ms), statistics.median(step_ms), max(step_ms)],
        "step_spread_50": ({"ms_min_p10_median_p90_max": [spread_ms[0], spread_ms[len(spread_ms) // 10],
                                                           statistics.median(spread_ms),
                                                           spread_ms[(9 * len(spread_ms)) // 10], spread_ms[-1]],
                            "us_per_layer_median": statistics.median(spread_ms) * 1e3 / st.L,
                            "note": "50 more graph replays after the timed region, each with its own queries"}
                           if spread_ms else None),
        "e2e_step_ms_min_median_max": [min(e2e_steps) * 1e3, statistics.median(e2e_steps) * 1e3,
                                       max(e2e_steps) * 1e3],
        "wall_ms_per_step": (wall1 - wall0) * 1e3 / args.steps,
        "eager_issue_us_per_layer": issue_s * 1e6 / st.L,
        "clocks": clk,
    }
    if hbm_scan is not None:
        line["hbm_scan"] = hbm_scan
    if fixed136 is not None:
        if "us_per_layer" in fixed136:
            fixed136["speedup_of_fathom"] = fixed136["us_per_layer"] / us_layer
            fixed136["note"] = ("the 32 channels of largest g at depth 4 (128 code bits + 8 scale bits per token) "
                                "through the same kernels and path; the pages report 1.67x at 1M tokens on an "
                                "A100 with PCIe 4.0 (Tab. 2), context only")
        line["vs_136bit"] = fixed136
    if st.host:
        line["link_gbs_peak"] = link_gbs
        line["link_gbs_sm_loads"] = sm_link_gbs
        line["link_roofline_frac_of_step"] = (scanned / (link_gbs * 1e9)) / (elapsed / (args.steps * L))
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.budget)
        try:
            line["cpu_baseline"]["all_cores"] = cpu_baseline_parallel(w, args.budget)
        except Exception as exc:   # reported as missing, never as a number
            log(f"[bench] all-cores CPU baseline unavailable: {exc}")
            line["cpu_baseline"]["all_cores"] = {"error": str(exc)[:200]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
