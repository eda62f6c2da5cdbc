"""The C-ABI library loads and exports every symbol include/fathom.h declares,
and argument validation rejects bad calls before any CUDA work (no GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

from bit_plane_kv_gb300 import binding as B
from bit_plane_kv_gb300 import build as BUILD

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fathom.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fathom_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    BUILD.build()
    return B.lib()


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert len(syms) >= 10, syms
    for s in syms:
        assert hasattr(lib, s), s
    # and the binding knows every one of them
    assert sorted(B.SIGNATURES) == syms


def test_version_and_struct_sizes(lib):
    assert "sm_103a" in B.version()
    assert ctypes.sizeof(B.Shape) == 9 * 4
    assert B.RUN_BYTES == 24


def rc_msg(lib, rc):
    return rc, lib.fathom_last_error().decode()


@pytest.mark.parametrize("field,value,frag", [
    ("units", 0, "units"), ("n", 0, "n must"), ("D", 0, "D must"), ("D", 129, "D must"),
    ("G", 3, "G must"), ("k", 0, "k must"), ("k", 5000, "k must"), ("n_sink", -1, "n_sink"),
    ("n_cap", 100, "n_cap"), ("scan_ctas_per_sm", -1, "scan_ctas_per_sm"), ("scan_ctas_per_sm", 9, "scan_ctas_per_sm"),
])
def test_shape_validation(lib, field, value, frag):
    s = B.make_shape(2, 4096, 128, 4, 64)
    setattr(s, field, value)
    dummy = ctypes.c_void_p(16)   # never dereferenced: validation fails first
    rc = lib.fathom_scan_topk(ctypes.byref(s), dummy, dummy, 0, 0, 0, dummy, dummy, dummy, dummy,
                              None, dummy, 1 << 30, None)
    rc, msg = rc_msg(lib, rc)
    assert rc == 1 and frag in msg, msg


def test_forced_exceeds_k(lib):
    s = B.make_shape(1, 4096, 128, 4, 20, 4, 32)
    assert lib.fathom_workspace_size(ctypes.byref(s), 0) == 0
    assert "forced" in lib.fathom_last_error().decode()


def test_null_pointers_and_small_workspace(lib):
    s = B.make_shape(1, 4096, 128, 4, 64)
    dummy = ctypes.c_void_p(256)
    rc = lib.fathom_quantize_pack(ctypes.byref(s), None, 0, dummy, dummy, None)
    assert rc_msg(lib, rc) == (1, "keys is NULL")
    need = lib.fathom_workspace_size(ctypes.byref(s), B.WS_SCAN_TOPK)
    assert need > 0
    rc = lib.fathom_scan_topk(ctypes.byref(s), dummy, dummy, 0, 0, 0, dummy, dummy, dummy, dummy,
                              None, dummy, need - 1, None)
    rc, msg = rc_msg(lib, rc)
    assert rc == 3 and "workspace too small" in msg
    rc = lib.fathom_scan_topk(ctypes.byref(s), dummy, dummy, 7, 0, 0, dummy, dummy, dummy, dummy,
                              None, dummy, need, None)
    assert rc_msg(lib, rc)[0] == 1
    rc = lib.fathom_plan_fixed(ctypes.byref(s), dummy, dummy, 0, 4, dummy, dummy, None)
    assert rc_msg(lib, rc)[0] == 1
    rc = lib.fathom_calibrate(1, 1, 128, dummy, None, dummy, None)
    assert rc_msg(lib, rc)[0] == 1
    rc = lib.fathom_sparse_attn(ctypes.byref(s), dummy, dummy, dummy, dummy, dummy, dummy,
                                lib.fathom_workspace_size(ctypes.byref(s), 1) - 1, None)
    assert rc_msg(lib, rc)[0] == 3


def test_workspace_sizes_scale_with_shape(lib):
    small = B.make_shape(1, 4096, 128, 4, 64)
    big = B.make_shape(8, 1 << 20, 128, 4, 512)
    assert 0 < B.workspace_size(small, 0) < B.workspace_size(big, 0)
    assert 0 < B.workspace_size(small, 1) <= B.workspace_size(big, 1)
    assert 0 < B.workspace_size(small, 2) <= B.workspace_size(big, 2)
    assert 0 < B.workspace_size(small, 3) <= B.workspace_size(big, 3)
    assert B.workspace_size(big, 4) == 0


def _attn_rows(pairs, k, sms=152):
    # kept-list entries per attention CTA for `pairs` grid rows of one head (the
    # library's rule; without a device it assumes 152 SMs)
    ctas128 = pairs * -(-k // 128)
    ctas512 = pairs * -(-k // 512)
    return 512 if ctas512 >= 4 * sms else (256 if ctas128 > 4 * sms else 128)


@pytest.mark.parametrize("units,G,k,D", [(1, 4, 64, 128), (8, 4, 512, 128), (39, 4, 512, 128), (152, 4, 512, 128),
                                         (256, 4, 512, 128), (16387, 4, 40, 128), (3, 8, 2048, 98), (5, 2, 300, 64)])
def test_attention_workspace_covers_both_launch_forms(lib, units, G, k, D):
    # the union form (one grid row per unit, G heads) and the per-head form (one grid
    # row per unit and head) share one workspace: partial states of whichever needs
    # more, then a ticket per (unit, head)
    shape = B.make_shape(units, 4096, D, G, k)
    ru = _attn_rows(units * G, k)                  # union form: units rows of G heads each
    rh = _attn_rows(units * G, k)                  # per-head form: units x G rows of one head
    splits_union = G * -(-k // ru)
    splits_head = -(-k // rh)
    part = max(units * splits_union * G, units * G * splits_head) * (D + 2) * 4
    align = lambda x: (x + 255) // 256 * 256
    need = align(align(part) + units * G * 4)
    assert B.workspace_size(shape, 1) == need


def test_fidelity_reference_calls_validate_arguments(lib):
    d = ctypes.c_void_p(256)
    s = B.make_shape(2, 4096, 128, 4, 64)
    need = lib.fathom_workspace_size(ctypes.byref(s), B.WS_SCAN_TOPK)
    rc = lib.fathom_exact_topk(ctypes.byref(s), None, d, d, d, None, d, need, None)
    assert rc_msg(lib, rc)[0] == 1
    rc = lib.fathom_exact_topk(ctypes.byref(s), d, d, d, d, None, d, need - 1, None)
    assert rc_msg(lib, rc)[0] == 3
    dn = lib.fathom_workspace_size(ctypes.byref(s), B.WS_DENSE_ATTN)
    rc = lib.fathom_dense_attn(ctypes.byref(s), d, d, d, None, d, dn, None)
    assert rc_msg(lib, rc) == (1, "out is NULL")
    rc = lib.fathom_dense_attn(ctypes.byref(s), d, d, d, d, d, dn - 1, None)
    assert rc_msg(lib, rc)[0] == 3


def test_rotated_basis_calls_validate_arguments(lib):
    d = ctypes.c_void_p(256)
    rc = lib.fathom_calibrate_klt(1, 1, 128, d, d, d, d, None)
    assert rc_msg(lib, rc)[0] == 1 and "m >= 2" in lib.fathom_last_error().decode()
    rc = lib.fathom_calibrate_klt(1, 16, 128, d, None, d, d, None)
    assert rc_msg(lib, rc) == (1, "mean is NULL")
    s = B.make_shape(2, 4096, 128, 4, 64)
    rc = lib.fathom_rotate_keys(ctypes.byref(s), d, 0, 0, d, d, d, None)
    assert rc_msg(lib, rc)[0] == 1 and "groups" in lib.fathom_last_error().decode()
    rc = lib.fathom_rotate_keys(ctypes.byref(s), d, 7, 1, d, d, d, None)
    assert rc_msg(lib, rc)[0] == 1
    rc = lib.fathom_rotate_query(ctypes.byref(s), d, 1, d, None, None)
    assert rc_msg(lib, rc) == (1, "q_rot is NULL")


def test_append_block_validates_its_block(lib):
    d = ctypes.c_void_p(256)
    s = B.make_shape(2, 4096, 128, 4, 64, n_cap=4160)
    for block, count in ((-1, 64), (0, 0), (0, 65), (65, 1), (64, 65)):
        rc = lib.fathom_append_block(ctypes.byref(s), d, 1, block, count, d, d, None)
        assert rc_msg(lib, rc)[0] == 1 and "append_block" in lib.fathom_last_error().decode()
    rc = lib.fathom_append_block(ctypes.byref(s), d, 1, 65, 0, d, d, None)
    assert rc_msg(lib, rc)[0] == 1


def test_online_basis_validates_arguments(lib):
    d = ctypes.c_void_p(256)
    s = B.make_shape(2, 4096, 128, 4, 64)
    need = lib.fathom_workspace_size(ctypes.byref(s), B.WS_KLT_ONLINE)
    assert need > 0
    rc = lib.fathom_klt_online(ctypes.byref(s), d, None, d, d, d, need, None)
    assert rc_msg(lib, rc) == (1, "mean is NULL")
    rc = lib.fathom_klt_online(ctypes.byref(s), d, d, d, d, d, need - 1, None)
    assert rc_msg(lib, rc)[0] == 3
    one = B.make_shape(2, 1, 128, 4, 1, 0, 0)
    rc = lib.fathom_klt_online(ctypes.byref(one), d, d, d, d, d, need, None)
    assert rc_msg(lib, rc)[0] == 1 and "n >= 2" in lib.fathom_last_error().decode()


def test_plane_key_attention_validates_arguments(lib):
    d = ctypes.c_void_p(256)
    s = B.make_shape(2, 4096, 128, 4, 64)
    need = lib.fathom_workspace_size(ctypes.byref(s), B.WS_SPARSE_ATTN)
    rc = lib.fathom_sparse_attn_planes(ctypes.byref(s), None, d, d, d, d, d, d, need, None)
    assert rc_msg(lib, rc) == (1, "planes is NULL")
    rc = lib.fathom_sparse_attn_planes(ctypes.byref(s), d, d, d, d, d, d, d, need - 1, None)
    assert rc_msg(lib, rc)[0] == 3


def test_fidelity_helpers_validate_and_greedy_matches_oracle(lib):
    # rows == 0 enqueues nothing; bad sizes are rejected before any launch
    assert lib.fathom_rel_err(0, 128, None, None, None, None) == 0
    assert rc_msg(lib, lib.fathom_rel_err(4, 0, None, None, None, None))[0] == 1
    assert rc_msg(lib, lib.fathom_set_overlap(4, 0, None, None, None, None))[0] == 1
    assert lib.fathom_set_overlap(0, 8, None, None, None, None) == 0
    # the greedy allocation is host code: it runs here and must equal the oracle's
    from oracle import oracle as O
    rng = np.random.default_rng(41)
    for trial in range(40):
        L, levels = int(rng.integers(1, 9)), int(rng.integers(1, 15))
        err = rng.uniform(0, 1, size=(L, levels))
        if trial % 3 == 0:
            err = np.round(err, 1)                        # many ties
        for b_mean in sorted({24, 24 + 8 * (levels - 1), 24 + 8 * int(rng.integers(0, levels))}):
            np.testing.assert_array_equal(B.fathom_greedy_budgets(err, 24, 8, b_mean),
                                          O.greedy_budgets(err, 24, 8, b_mean))
    with pytest.raises(B.FathomError):
        B.fathom_greedy_budgets(np.zeros((2, 14)), 24, 8, 50)           # 50 is not a level
    with pytest.raises(B.FathomError):
        B.fathom_greedy_budgets(np.full((2, 14), np.nan), 24, 8, 48)
    with pytest.raises(B.FathomError):
        B.fathom_greedy_budgets(np.zeros((2, 3)), 24, 8, 48)            # above the top level (40)


def test_debug_status_reports_a_build_without_checks(lib):
    # the default build compiles every bounds check away: the call says so and writes zeros
    out = (ctypes.c_uint64 * 3)(7, 7, 7)
    rc = lib.fathom_debug_status(0, ctypes.cast(out, ctypes.c_void_p))
    code, msg = rc_msg(lib, rc)
    assert code == 1 and "without the debug checks" in msg
    assert list(out) == [0, 0, 0]
    assert rc_msg(lib, lib.fathom_debug_status(3, ctypes.cast(out, ctypes.c_void_p)))[0] == 1
    assert rc_msg(lib, lib.fathom_debug_status(0, None)) == (1, "first_failure is NULL")


# ---- the scan's grid choice, seen through the workspace size (host logic, no device:
# the library then assumes 152 SMs with 3 resident scan CTAs each)
def _scan_makespan(units, n_sub, chunks, slots, unit_fast):
    import heapq
    total = units * chunks
    ctr = [0] * units
    took = [False] * total
    q = [(0.0, i) for i in range(min(total, slots))]
    heapq.heapify(q)
    nxt, end = min(total, slots), 0.0
    while q:
        t, i = heapq.heappop(q)
        u = i % units if unit_fast else i // chunks
        if ctr[u] < n_sub:
            ctr[u] += 1
            took[i] = True
            heapq.heappush(q, (t + 1.0, i))
            continue
        t2 = t + (1.0 if took[i] else 0.1)
        end = max(end, t2)
        if nxt < total:
            heapq.heappush(q, (t2, nxt))
            nxt += 1
    return end


def _scan_chunks(units, n, slots=152 * 3):
    n_sub = -(-(-(-n // 64)) // 32)
    best, best_cost = 1, None
    for c in range(1, min(n_sub, 4096) + 1):
        waves = -(-(units * c) // slots)
        cost = waves * (-(-n_sub // c) + 1)
        if best_cost is None or cost < best_cost:
            best, best_cost = c, cost
        if units * c >= 8 * slots:
            break
    if units < slots and slots % units and units * n_sub <= 1000000:
        q0 = slots // units + 1
        uf_cost, uf_best = best_cost, 0
        for c in range(q0, min(4 * q0, n_sub, 4096) + 1):
            t = _scan_makespan(units, n_sub, c, slots, True)
            if t < uf_cost:
                uf_cost, uf_best = t, c
        if uf_best:
            best = uf_best
    return best


def _scan_ws(units, n, G, k, chunks, n_sink=4, n_recent=32):
    a = lambda x: (x + 255) // 256 * 256
    ns = min(n_sink, n)
    r0 = max(ns, n - n_recent)
    nf = ns + n - r0
    ksel = max(k - nf, 0)
    cap = a(ksel + 256 + 2 * 2048)
    ks1 = max(ksel, 1)
    m = min(max(-(-4 * ks1 // chunks), 32), ks1)
    parts = max(min(-(-(chunks * 3 * m) // 8192), chunks, 1024), 1)
    ctas, uh = units * chunks, units * G
    off = a(ctas * G * cap * 8)
    off = a(off + ctas * G * 4)
    off = a(off + ctas * G * 8)
    off = a(off + ctas * G * 4)
    off = a(off + uh * max(nf, 1) * 4)
    off = a(off + uh * parts * ks1 * 8)
    off = a(off + uh * parts * 4)
    off = a(off + uh * 4)
    off = a(off + uh * 4)
    n_sub = -(-(-(-n // 64)) // 32)
    off = a(off + units * 4)
    return a(off + units * n_sub * 4)


@pytest.mark.parametrize("units,n", [(8, 1 << 20), (8, 1 << 15), (256, 1 << 16), (300, 1 << 16), (100, 1 << 17),
                                     (2048, 1 << 16), (1, 4096), (24, 1 << 20)])
def test_scan_grid_choice_matches_a_simulation_of_the_schedule(lib, units, n):
    # the chunk count behind the workspace size is the one a direct simulation of
    # the shared sub-chunk counters picks (unit-fastest launch only where the units
    # do not fill the resident slots evenly); for 256 units of 64k tokens it is the
    # unit-fastest launch with 8 CTAs per unit
    G, k = 4, 512
    shape = B.make_shape(units, n, 128, G, k)
    got = B.workspace_size(shape, 0)
    c = _scan_chunks(units, n)
    assert got == _scan_ws(units, n, G, k, c), (units, n, c)
    if (units, n) == (256, 1 << 16):
        assert c == 8
